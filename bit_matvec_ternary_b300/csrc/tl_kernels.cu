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
//   Work.  The launch's (16-row tile, 128-column block) units are ordered row
//   tile by row tile; CTA c owns the contiguous range [c*Lc, (c+1)*Lc), so
//   every CTA streams the same number of bytes and a row tile spans at most
//   two CTAs.  Inside a CTA the k-range is processed in passes of KS blocks
//   (the activations of one pass fit the staging buffer at 8 tokens); the 16
//   warps split each pass's units into contiguous ranges.
//   Weights.  Each warp streams its units with cp.async.bulk into its own
//   ring of shared-memory slots (up to 4 tiles, 2 KB, per copy, completing
//   on the slot's mbarrier), running ahead across passes.  A TL2P v1 tile is
//   in mma.m16n8k16 A-fragment order: register f of a 16-column step is
//   (word << 2q) & 0xC000C000, a bf16x2 pair of +-2.0 / +-0.0 -- one shift
//   (IMAD, FMA pipe) and one AND (LOP3, ALU pipe) per two weights; the
//   tensor cores do the multiply-adds (products exact, fp32 sums).
//   Activations.  Staged per pass in shared memory in B-fragment order (mode
//   B converts int8 to bf16, exact); columns n >= N repeat token N-1 and
//   their results are discarded, so no lane is predicated off.
//   Reduction.  A warp that covers all of a row tile's units in a pass adds
//   its sum straight into the CTA's row accumulator (shared memory); rows
//   split between warps go through per-warp boundary slots that are added in
//   warp order after the pass.  A row tile cut by a CTA boundary is finished
//   by whichever of its two CTAs arrives second (workspace counter), adding
//   the two halves in a fixed order.  The plan never depends on N, so every
//   token's result is bitwise independent of the batch.

#include "tl.h"
#include "tl_internal.cuh"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <algorithm>
#include <cstring>

namespace {

constexpr int kWarps = 16;            // warps per CTA of the N <= 8 kernel (one CTA per SM)
constexpr int kThreads = kWarps * 32;
constexpr int kChunkTiles = 4;        // tiles (512 B each) per bulk copy
constexpr int kSlots = 2;             // bulk copies in flight per warp
constexpr int kRingBytes = kWarps * kSlots * kChunkTiles * 512;   // 64 KB
constexpr int kNMax = 8;              // tokens per launch (mma n = 8)
constexpr int kMaxDevices = 64;
constexpr int kStageBlocks = 16;      // 128-column blocks per pass (32 KB at 8 tokens)
constexpr int kMaxCtaRows = 32;       // row tiles one CTA may touch
constexpr long long kWaitLimit = 1ll << 31;   // SM cycles before a wait gives up

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
    int KS;         // blocks per pass
    int S;          // passes
    int K;
    int U;          // units = R * KB
    int Lc;         // units per CTA (the last CTAs may get fewer)
    const void *X;  // bf16 [N][K] (mode A) or int8 [N][K] (mode B)
    const float *s;
    const int32_t *z;
    int N;
    int mode;
    int out;
    float *part;    // halves of CTA-split row tiles [R][2][N][16]
    unsigned long long *cnt;  // [R] blocks arrived; zero between launches
    int *status;    // workspace status word
};

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
// The CTA's unit range and the row tiles it touches.
struct CtaGeo {
    int cu0, cu1;           // units [cu0, cu1), unit = row_tile * KB + block
    int r_first, r_last;    // row tiles touched (r_last < r_first: none)
    int lo_first, hi_last;  // first block of r_first, one past the last block of r_last
};

__device__ __forceinline__ CtaGeo cta_geo(const GroupArgs &a, int c) {
    CtaGeo g;
    g.cu0 = min(c * a.Lc, a.U);
    g.cu1 = min(g.cu0 + a.Lc, a.U);
    if (g.cu1 > g.cu0) {
        g.r_first = g.cu0 / a.KB;
        g.r_last = (g.cu1 - 1) / a.KB;
        g.lo_first = g.cu0 - g.r_first * a.KB;
        g.hi_last = g.cu1 - g.r_last * a.KB;
    } else {
        g.r_first = 0; g.r_last = -1; g.lo_first = 0; g.hi_last = 0;
    }
    return g;
}

// Blocks [lo, hi) of row tile r that the CTA covers in pass s.
__device__ __forceinline__ void row_span(const GroupArgs &a, const CtaGeo &g, int r, int s,
                                         int &lo, int &hi) {
    lo = max(r == g.r_first ? g.lo_first : 0, s * a.KS);
    hi = min(r == g.r_last ? g.hi_last : a.KB, (s + 1) * a.KS);
}

__device__ __forceinline__ int row_count(const GroupArgs &a, const CtaGeo &g, int r, int s) {
    int lo, hi;
    row_span(a, g, r, s, lo, hi);
    return max(0, hi - lo);
}

__device__ __forceinline__ int pass_units(const GroupArgs &a, const CtaGeo &g, int s) {
    if (g.r_last < g.r_first) return 0;
    const int c0 = row_count(a, g, g.r_first, s);
    if (g.r_last == g.r_first) return c0;
    return c0 + (g.r_last - g.r_first - 1) * a.KS + row_count(a, g, g.r_last, s);
}

// Row tile and block of the i-th unit of pass s in the CTA.
__device__ __forceinline__ void pass_locate(const GroupArgs &a, const CtaGeo &g, int s, int i,
                                            int &r, int &b) {
    int lo, hi;
    row_span(a, g, g.r_first, s, lo, hi);
    const int c0 = max(0, hi - lo);
    if (i < c0) { r = g.r_first; b = lo + i; return; }
    const int j = i - c0;
    const int mid = g.r_last > g.r_first ? (g.r_last - g.r_first - 1) * a.KS : 0;
    if (j < mid) { r = g.r_first + 1 + j / a.KS; b = s * a.KS + j % a.KS; return; }
    row_span(a, g, g.r_last, s, lo, hi);
    r = g.r_last;
    b = lo + (j - mid);
}

// A warp's walk over its units, pass after pass, in chunks: runs of at most
// kChunkTiles consecutive blocks of one row tile (contiguous in memory).
struct Walk {
    int s, i, iend;          // pass, unit index in the pass, end of the warp's range
    int r, b, row_hi;        // current row tile, block, end block of the row in this pass
    int gi, rl;              // matrix of the group and its local row tile
    int n;                   // tiles in the current chunk (0: done)

    __device__ void map_row(const GroupArgs &a) {
        gi = 0;
        while (gi + 1 < a.G && a.rt_off[gi + 1] <= r) ++gi;
        rl = r - a.rt_off[gi];
    }
    __device__ void enter(const GroupArgs &a, const CtaGeo &g, int w) {
        // from pass s on: the first pass in which warp w has units
        for (; s < a.S; ++s) {
            const int np = pass_units(a, g, s);
            const int lw = (np + kWarps - 1) / kWarps;
            i = min(w * lw, np);
            iend = min(i + lw, np);
            if (i < iend) {
                pass_locate(a, g, s, i, r, b);
                int lo;
                row_span(a, g, r, s, lo, row_hi);
                map_row(a);
                n = min(kChunkTiles, min(iend - i, row_hi - b));
                return;
            }
        }
        n = 0;
    }
    __device__ void start(const GroupArgs &a, const CtaGeo &g, int w) {
        s = 0;
        enter(a, g, w);
    }
    __device__ void next(const GroupArgs &a, const CtaGeo &g, int w) {
        i += n;
        b += n;
        if (i >= iend) {
            ++s;
            enter(a, g, w);
            return;
        }
        if (b >= row_hi) {
            ++r;
            int lo;
            row_span(a, g, r, s, lo, row_hi);
            b = lo;
            map_row(a);
        }
        n = min(kChunkTiles, min(iend - i, row_hi - b));
    }
    __device__ __forceinline__ const char *src(const GroupArgs &a) const {
        return a.packed[gi] + ((long long)rl * a.KB + b) * 512;
    }
};

// ------------------------------------------------------------ epilogue
// Y[n][m] from acc_y = sum_k w*x (mode A) or the exact integer sum_k w*q (mode B).
__device__ __forceinline__ void store_out(const GroupArgs &a, int gi, int m, int n, float acc) {
    const int M = a.M[gi];
    float y;
    if (a.mode == TL_MODE_BF16) {
        y = __fmul_rn(acc, a.scale[gi][m]);
    } else {
        const int iacc = __float2int_rn(acc);
        if (a.out == TL_OUT_I32_RAW) {
            reinterpret_cast<int32_t *>(a.Y[gi])[(long long)n * M + m] = iacc;
            return;
        }
        const int corrected = iacc - a.z[n] * a.rowsum[gi][m];
        y = __fmul_rn(__fmul_rn((float)corrected, a.s[n]), a.scale[gi][m]);
    }
    if (a.out == TL_OUT_F32)
        reinterpret_cast<float *>(a.Y[gi])[(long long)n * M + m] = y;
    else
        reinterpret_cast<__nv_bfloat16 *>(a.Y[gi])[(long long)n * M + m] = __float2bfloat16_rn(y);
}

// The 16 x N results of row tile r held as acc[n * 16 + row] (sums of +-2
// weights: halved here, exactly).  One warp; lane (g, t) stores rows g, g+8
// of tokens 2t, 2t+1.
__device__ __forceinline__ void store_row_tile(const GroupArgs &a, int r, const float *acc,
                                               int lane) {
    const int g = lane >> 2, t = lane & 3;
    int gi = 0;
    while (gi + 1 < a.G && a.rt_off[gi + 1] <= r) ++gi;
    const int rl = r - a.rt_off[gi];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int m = rl * 16 + g + 8 * h, n = 2 * t + e;
            if (m < a.M[gi] && n < a.N) store_out(a, gi, m, n, acc[n * 16 + g + 8 * h] * 0.5f);
        }
}

// One 128-column block of one 16-row tile: 8 MMAs over the lane's 16-byte
// slice of the tile (w) and the 4 B-fragment quarters (b).
__device__ __forceinline__ void tile_mma(float (&c)[4][4], const uint4 &w, const uint4 (&b)[4]) {
    const uint32_t M2 = 0xC000C000u;
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
    // four independent accumulator chains; consecutive MMAs never share one
#pragma unroll
    for (int qd = 0; qd < 4; ++qd)
        mma_bf16_16816(c[qd], wd[qd] & M2, (wd[qd] << 2) & M2, (wd[qd] << 4) & M2,
                       (wd[qd] << 6) & M2, b[qd].x, b[qd].y);
#pragma unroll
    for (int qd = 0; qd < 4; ++qd)
        mma_bf16_16816(c[qd], (wd[qd] << 8) & M2, (wd[qd] << 10) & M2, (wd[qd] << 12) & M2,
                       (wd[qd] << 14) & M2, b[qd].z, b[qd].w);
}

// ------------------------------------------------------------ kernel
// kModeA: bf16 activations (else int8 from the quantiser).  NT: token
// columns staged (a power of two >= N).
template <bool kModeA, int NT>
__global__ void __launch_bounds__(kThreads)
tl_mma_kernel(const __grid_constant__ GroupArgs a) {
    constexpr int XQ = NT * 4;                  // uint4 per 32-column quarter
    constexpr int XB = 4 * XQ;                  // uint4 per 128-column block
    constexpr int RV = 16 * NT;                 // floats per row-tile result
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;                                              // [kWarps][kSlots][2 KB]
    uint4 *xs = reinterpret_cast<uint4 *>(smem + kRingBytes);          // one pass of X
    float *acc = reinterpret_cast<float *>(smem + kRingBytes + a.KS * XB * 16);  // [rows][RV]
    __shared__ float bslot[kWarps][2][RV];      // boundary pieces of the current pass
    __shared__ int bslot_row[kWarps][2];
    __shared__ __align__(8) unsigned long long bars[kWarps][kSlots];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const CtaGeo geo = cta_geo(a, blockIdx.x);
    const int nrows = geo.r_last - geo.r_first + 1;
    const int N = a.N;

    if (threadIdx.x < kWarps * kSlots)
        mbar_init(smem_u32(&bars[0][0]) + 8u * threadIdx.x, 1);
    if (threadIdx.x < kWarps * 2) (&bslot_row[0][0])[threadIdx.x] = -1;
    for (int i = threadIdx.x; i < nrows * RV; i += kThreads) acc[i] = 0.f;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();

    // Weights do not depend on the previous kernel: start the bulk copies
    // before waiting for it.  The producer (lane 0) runs kSlots chunks ahead
    // of the consumer, across pass boundaries.
    const uint32_t ring_w = smem_u32(ring) + warp * (kSlots * kChunkTiles * 512);
    const uint32_t bar_w = smem_u32(&bars[warp][0]);
    Walk pf;
    pf.start(a, geo, warp);
    if (lane == 0)
        for (int k = 0; k < kSlots && pf.n > 0; ++k) {
            bulk_load(ring_w + k * (kChunkTiles * 512), pf.src(a), pf.n * 512, bar_w + 8u * k);
            pf.next(a, geo, warp);
        }
    griddep_wait();
    griddep_launch();

    Walk cw;
    cw.start(a, geo, warp);
    int slot = 0;
    uint32_t phases = 0;                        // parity bit per slot
    bool ok = true;
    float c[4][4];

    for (int s = 0; s < a.S; ++s) {
        // ---- stage X for pass s in B-fragment order:
        // word ((((bp*4 + qd)*NT + n)*4 + t)*4 + w) holds x[n'][k], x[n'][k+1],
        // n' = min(n, N-1), k = (s*KS + bp)*128 + 16*(2qd + w/2) + 2t + 8*(w%2).
        {
            const int words = a.KS * 64 * NT;
            uint32_t *xw = reinterpret_cast<uint32_t *>(xs);
            for (int idx = threadIdx.x; idx < words; idx += kThreads) {
                const int w = idx & 3, tt = (idx >> 2) & 3;
                const int n = min((idx >> 4) % NT, N - 1);
                const int rest = (idx >> 4) / NT;
                const int qd = rest & 3, bp = rest >> 2;
                const int k = (s * a.KS + bp) * 128 + 16 * (2 * qd + (w >> 1)) + 2 * tt + 8 * (w & 1);
                uint32_t lo = 0, hi = 0;
                if (kModeA) {
                    const uint16_t *x = reinterpret_cast<const uint16_t *>(a.X) + (long long)n * a.K;
                    if (k < a.K) lo = x[k];
                    if (k + 1 < a.K) hi = x[k + 1];
                } else {
                    const int8_t *x = reinterpret_cast<const int8_t *>(a.X) + (long long)n * a.K;
                    if (k < a.K) lo = __bfloat16_as_ushort(__float2bfloat16_rn((float)x[k]));
                    if (k + 1 < a.K) hi = __bfloat16_as_ushort(__float2bfloat16_rn((float)x[k + 1]));
                }
                xw[idx] = lo | (hi << 16);
            }
        }
        __syncthreads();

        // ---- this warp's units of pass s
        int run_lo = cw.b, nslot = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
        while (ok && cw.n > 0 && cw.s == s) {
            const bool got = __all_sync(0xffffffffu,
                                        mbar_wait(bar_w + 8u * slot, (phases >> slot) & 1u, a.status));
            if (!got) { ok = false; break; }
            phases ^= 1u << slot;
            const uint4 *tiles = reinterpret_cast<const uint4 *>(
                ring + warp * (kSlots * kChunkTiles * 512) + slot * (kChunkTiles * 512)) + lane;
            const uint4 *xb = xs + (cw.b - s * a.KS) * XB + (g % NT) * 4 + t;
            if (cw.n == kChunkTiles) {
                // full chunk: load tile i+1 while tile i is multiplied
                uint4 w = tiles[0];
                uint4 bq[4];
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) bq[qd] = xb[qd * XQ];
#pragma unroll
                for (int i = 0; i < kChunkTiles; ++i) {
                    uint4 wn = w, bn[4] = {bq[0], bq[1], bq[2], bq[3]};
                    if (i + 1 < kChunkTiles) {
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
                for (int i = 0; i < cw.n; ++i) {
                    const uint4 w = tiles[i * 32];
                    uint4 bq[4];
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd) bq[qd] = xb[i * XB + qd * XQ];
                    tile_mma(c, w, bq);
                }
            }
            // end of a run of one row tile: this chunk ends the row or the warp's range
            const bool run_end = (cw.b + cw.n == cw.row_hi) || (cw.i + cw.n == cw.iend);
            if (run_end) {
                float v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) v[q] = (c[0][q] + c[1][q]) + (c[2][q] + c[3][q]);
                int lo, hi;
                row_span(a, geo, cw.r, s, lo, hi);
                const int rho = cw.r - geo.r_first;
                // lane (g, t) holds rows g, g+8 of tokens 2t, 2t+1
                if (run_lo == lo && cw.b + cw.n == hi) {
                    // the whole row tile of this pass: no other warp touches it
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
                run_lo = cw.b + cw.n < cw.row_hi ? cw.b + cw.n : -1;   // next run starts a row
            }
            // refill this slot with the chunk kSlots ahead
            __syncwarp();
            if (lane == 0 && pf.n > 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                bulk_load(ring_w + slot * (kChunkTiles * 512), pf.src(a), pf.n * 512, bar_w + 8u * slot);
                pf.next(a, geo, warp);
            }
            cw.next(a, geo, warp);
            if (run_lo < 0) run_lo = cw.b;
            slot = slot + 1 == kSlots ? 0 : slot + 1;
        }
        __syncthreads();
        // ---- boundary pieces of pass s, added in warp order (one thread per element)
        if (threadIdx.x < RV) {
            for (int w = 0; w < kWarps; ++w)
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int rho = bslot_row[w][k];
                    if (rho >= 0) acc[rho * RV + threadIdx.x] += bslot[w][k][threadIdx.x];
                }
        }
        __syncthreads();
        if (threadIdx.x < kWarps * 2) (&bslot_row[0][0])[threadIdx.x] = -1;
        // (the next pass's staging __syncthreads orders this reset before reuse)
    }
    if (!ok) {
        // a copy never landed: drain what is still in flight (bounded), then leave
        for (int k = 0; k < kSlots; ++k) mbar_wait(bar_w + 8u * k, (phases >> k) & 1u, a.status);
        return;
    }

    // ---- results: rows covered entirely by this CTA go straight to Y; a row
    // tile cut by a CTA boundary is finished by the second of its two CTAs.
    for (int rho = warp; rho < nrows; rho += kWarps) {
        const int r = geo.r_first + rho;
        const int lo = r == geo.r_first ? geo.lo_first : 0;
        const int hi = r == geo.r_last ? geo.hi_last : a.KB;
        const float *v = acc + rho * RV;
        if (lo == 0 && hi == a.KB) {
            store_row_tile(a, r, v, lane);
            continue;
        }
        const int half = lo == 0 ? 0 : 1;       // 0: holds block 0 of the row
        float *dst = a.part + ((long long)r * 2 + half) * N * 16;
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
            const float *h0 = a.part + (long long)r * 2 * N * 16;
            // combine the halves (block-0 half first) through this CTA's acc row
            for (int e = lane; e < N * 16; e += 32)
                acc[rho * RV + e] = __ldcg(h0 + e) + __ldcg(h0 + N * 16 + e);
            __syncwarp();
            store_row_tile(a, r, acc + rho * RV, lane);
            if (lane == 0) a.cnt[r] = 0ull;
        }
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

constexpr int kMaxDynSmem = kRingBytes + kStageBlocks * 128 * kNMax * 2 + kMaxCtaRows * 16 * kNMax * 4;

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
                                             kMaxDynSmem) != cudaSuccess)
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
    int R, KB, KS, S, P, Lc, rows;
    long long U;
    size_t smem;       // dynamic shared memory for the given N
    size_t ws_bytes;   // workspace for the given N
};

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// The plan depends on the shapes and the SM count only, never on N, so every
// token is summed in the same order whatever the batch.
tl_status make_plan(const int *Ms, int G, int K, int N, int sms, Plan *p) {
    p->R = 0;
    for (int g = 0; g < G; ++g) p->R += (int)ceil_div(Ms[g], 16);
    p->KB = (int)ceil_div(K, 128);
    p->U = (long long)p->R * p->KB;
    if (p->U >= (1ll << 30)) return TL_ERR_SHAPE;
    // passes: the largest divisor of KB not above kStageBlocks
    p->KS = 1;
    for (int d = 1; d <= std::min(p->KB, kStageBlocks); ++d)
        if (p->KB % d == 0) p->KS = d;
    p->S = p->KB / p->KS;
    // CTAs: at most one per SM, and ranges of at least KB - 1 units so a row
    // tile never spans more than two CTAs
    long long P = sms;
    if (p->KB > 1) P = std::min<long long>(P, std::max<long long>(1, p->U / (p->KB - 1)));
    else P = std::min<long long>(P, p->U);
    p->P = (int)std::max<long long>(1, P);
    p->Lc = (int)ceil_div(p->U, p->P);
    p->rows = (int)(ceil_div(p->Lc + p->KB - 1, p->KB) + 1);
    p->rows = std::min(p->rows, p->R);
    if (p->rows > kMaxCtaRows) return TL_ERR_SHAPE;
    const int nt = padded_tokens(std::min(std::max(N, 1), kNMax));
    const int n = std::min(std::max(N, 1), kNMax);
    p->smem = (size_t)kRingBytes + (size_t)p->KS * 128 * nt * 2 + (size_t)p->rows * 16 * nt * 4;
    const size_t cnt_bytes = ((size_t)p->R * 8 + 255) / 256 * 256;
    p->ws_bytes = tl_internal::kStatusBytes + cnt_bytes + (size_t)p->R * 2 * 16 * n * 4;
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
        if (w.layout != TL_LAYOUT_TL2P_V1) return TL_ERR_UNSUPPORTED;
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
        return std::max(tl_internal::prefill_workspace_bytes(N, K, TL_MODE_BF16),
                        tl_internal::prefill_workspace_bytes(N, K, TL_MODE_I8));
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
    a.R = p.R; a.KB = p.KB; a.KS = p.KS; a.S = p.S; a.K = K; a.U = (int)p.U; a.Lc = p.Lc;
    const size_t xsz = mode == TL_MODE_BF16 ? 2 : 1;
    a.X = static_cast<const char *>(X) + (size_t)n0 * K * xsz;
    a.s = s ? s + n0 : nullptr;
    a.z = z ? z + n0 : nullptr;
    a.N = n; a.mode = mode; a.out = out;
    const size_t cnt_bytes = ((size_t)p.R * 8 + 255) / 256 * 256;
    char *wsb = static_cast<char *>(ws) + tl_internal::kStatusBytes;
    a.cnt = reinterpret_cast<unsigned long long *>(wsb);
    a.part = reinterpret_cast<float *>(wsb + cnt_bytes);
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
    *zeroed = kStatusBytes + ((size_t)p.R * 8 + 255) / 256 * 256;
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
