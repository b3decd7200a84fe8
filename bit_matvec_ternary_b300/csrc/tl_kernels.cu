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
//   Weights.  Each warp owns a contiguous range of (slice, 16-row tile,
//   128-column block) units and streams them with cp.async.bulk into its own
//   ring of shared-memory slots (one bulk copy moves up to 4 tiles, 2 KB,
//   and completes on the slot's mbarrier).  A TL2P v1 tile is in
//   mma.m16n8k16 A-fragment order: a lane's 16 bytes are 4 words, each
//   covering two 16-column steps, and register f of a step is
//   (word << 2q) & 0xC000C000, a bf16x2 pair of +-2.0 / +-0.0 -- one shift
//   (IMAD, FMA pipe) and one AND (LOP3, ALU pipe) per two weights.  The
//   tensor cores do the multiply-adds (bf16 x bf16 -> fp32, products exact).
//   Activations.  Staged once per CTA in shared memory in B-fragment order
//   (mode B converts int8 to bf16, exact).  Token columns n >= N read token
//   N-1 (their results are discarded), so no lane is predicated off.
//   Split-K.  Warp v owns units [v*L, min((v+1)*L, U)), L = ceil(U / warps).
//   A row tile whose k-range spans several warps is finished by the warp
//   that completes its arrival count (workspace counter); it adds the pieces
//   in a fixed order, so results are deterministic and every token's result
//   is independent of N.

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
constexpr int kSlots = 3;             // bulk copies in flight per warp
constexpr int kRingBytes = kWarps * kSlots * kChunkTiles * 512;   // 96 KB
constexpr int kNMax = 8;              // tokens per launch (mma n = 8)
constexpr int kMaxDevices = 64;
constexpr size_t kSmemLimit = 120 * 1024;   // activation staging budget per CTA
constexpr int kMaxSlice = 32;         // 128-column blocks per split-K slice, at most
constexpr int kMaxPending = 8;        // partial pieces a warp holds before publishing
constexpr int kMaxSlices = 32;        // split-K slices per launch (one flag bit each)
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
    int KS;         // blocks per slice
    int S;          // slices
    int K;
    long long U;    // units = R * KB
    long long V;    // warps in the grid
    int L;          // units per warp (the last warps may get fewer or none)
    const void *X;  // bf16 [N][K] (mode A) or int8 [N][K] (mode B)
    const float *s;
    const int32_t *z;
    int N;
    int mode;
    int out;
    float *part;    // split-K partials [R*S*2][N][16]
    unsigned long long *cnt;  // [R] arrivals: low 32 bits = blocks summed so far,
                              // bit 32+s = slice s arrived in two pieces; zero between launches
    int *status;    // workspace status word
};

__device__ __forceinline__ int bnd(const GroupArgs &a, int v) {
    return (int)min((long long)v * a.L, a.U);
}

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
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
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

// A run of consecutive tiles of one (slice, row tile) segment: at most
// kChunkTiles, never across a segment or the warp's range end, so its bytes
// are contiguous in the packed matrix.
struct Chunk {
    int u, s, r, bp, gi, rl, n;

    __device__ void seek(const GroupArgs &a, int u0, int u1) {
        u = u0;
        const int su = a.R * a.KS;
        s = u0 / su;
        const int rem = u0 - s * su;
        r = rem / a.KS;
        bp = rem - r * a.KS;
        gi = 0;
        while (gi + 1 < a.G && a.rt_off[gi + 1] <= r) ++gi;
        rl = r - a.rt_off[gi];
        size(a, u1);
    }
    __device__ __forceinline__ void size(const GroupArgs &a, int u1) {
        n = min(kChunkTiles, min(a.KS - bp, u1 - u));
    }
    __device__ __forceinline__ void next(const GroupArgs &a, int u1) {
        u += n;
        bp += n;
        if (bp == a.KS) {
            bp = 0;
            if (++r == a.R) {
                r = 0; ++s; gi = 0; rl = 0;
            } else if (r == a.rt_off[gi + 1]) {
                ++gi; rl = 0;
            } else {
                ++rl;
            }
        }
        size(a, u1);
    }
    __device__ __forceinline__ const char *src(const GroupArgs &a) const {
        return a.packed[gi] + ((long long)rl * a.KB + (long long)s * a.KS + bp) * 512;
    }
    __device__ __forceinline__ bool seg_end(const GroupArgs &a, int u1) const {
        return bp + n == a.KS || u + n == u1;
    }
};

// Y[n][m] from the scaled sum y_acc = sum_k w*x (mode A) or the exact
// integer sum_k w*q (mode B).
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

__device__ __forceinline__ void epilogue(const GroupArgs &a, int gi, int rl, int g, int t,
                                         const float (&c)[4]) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int m = rl * 16 + g + 8 * h;
            const int n = 2 * t + e;
            if (m < a.M[gi] && n < a.N) store_out(a, gi, m, n, c[2 * h + e]);
        }
}

// Sum every piece of row tile r in fixed (slice, piece) order and store Y.
// Called by the warp whose arrival completed the row tile's count; `split`
// has bit s set when slice s came in two pieces.
__device__ __noinline__ void reduce_row_tile(const GroupArgs &a, int r, unsigned split,
                                             int lane) {
    const int g = lane >> 2, t = lane & 3;
    int gi = 0;
    while (gi + 1 < a.G && a.rt_off[gi + 1] <= r) ++gi;
    const int rl = r - a.rt_off[gi];
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int ss = 0; ss < a.S; ++ss) {
        const int pieces = ((split >> ss) & 1u) ? 2 : 1;
        for (int pp = 0; pp < pieces; ++pp) {
            const float *src = a.part + (((long long)r * a.S + ss) * 2 + pp) * a.N * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int n = 2 * t + e;
                    if (n < a.N) acc[2 * h + e] += __ldcg(src + n * 16 + g + 8 * h);
                }
        }
    }
    epilogue(a, gi, rl, g, t, acc);
    if (lane == 0) a.cnt[r] = 0ull;
}

// Publish this warp's pending pieces.  The lanes' partial-sum stores are
// ordered before lane 0's counter update by __syncwarp, and the update is a
// release (and acquire) at GPU scope, so the warp that completes a row tile's
// count sees every piece; it then reduces the row tile.  No full fence.
__device__ __forceinline__ unsigned long long atomic_add_acq_rel(unsigned long long *p,
                                                                 unsigned long long v) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;"
                 : "=l"(old)
                 : "l"(p), "l"(v)
                 : "memory");
    return old;
}

__device__ __noinline__ void commit_pieces(const GroupArgs &a, const int *pend_r,
                                           const unsigned long long *pend_add, int count,
                                           int lane) {
    __syncwarp();
    for (int i = 0; i < count; ++i) {
        const int r = pend_r[i];
        unsigned long long now = 0ull;
        if (lane == 0) now = atomic_add_acq_rel(a.cnt + r, pend_add[i]) + pend_add[i];
        now = __shfl_sync(0xffffffffu, now, 0);
        if ((unsigned)(now & 0xffffffffull) == (unsigned)a.KB) {
            __syncwarp();
            reduce_row_tile(a, r, (unsigned)(now >> 32), lane);
        }
    }
}

// Emit one piece (row tile r, slice s, piece p, nk blocks): the final result
// when it covers the whole k-range, else its partial sums go to the workspace
// and the piece joins the warp's pending list.  Returns the new list length.
__device__ __noinline__ int emit_piece(const GroupArgs &a, int r, int s, int p, int nk, int gi,
                                       int rl, int lane, float c0, float c1, float c2, float c3,
                                       int *pend_r, unsigned long long *pend_add,
                                       int pend_count) {
    const int g = lane >> 2, t = lane & 3;
    const float c[4] = {c0, c1, c2, c3};
    if (a.S == 1 && nk == a.KB) {   // the whole k-range in one piece: final
        epilogue(a, gi, rl, g, t, c);
        return pend_count;
    }
    const long long slot = ((long long)r * a.S + s) * 2 + p;
    float *dst = a.part + slot * a.N * 16;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = 2 * t + e;
            if (n < a.N) __stcg(dst + n * 16 + g + 8 * h, c[2 * h + e]);
        }
    if (lane == 0) {
        pend_r[pend_count] = r;
        pend_add[pend_count] = (unsigned long long)nk | ((unsigned long long)p << (32 + s));
    }
    __syncwarp();
    if (++pend_count == kMaxPending) {
        commit_pieces(a, pend_r, pend_add, pend_count, lane);
        pend_count = 0;
    }
    return pend_count;
}

// One 128-column block of one 16-row tile: 8 MMAs over the lane's 16-byte
// slice of the tile (w) and the 4 B-fragment quarters (b).
__device__ __forceinline__ void tile_mma(float (&c)[4][4], const uint4 &w, const uint4 (&b)[4]) {
    const uint32_t M2 = 0xC000C000u;
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
        const uint32_t word = qd == 0 ? w.x : qd == 1 ? w.y : qd == 2 ? w.z : w.w;
        mma_bf16_16816(c[qd], word & M2, (word << 2) & M2, (word << 4) & M2, (word << 6) & M2,
                       b[qd].x, b[qd].y);
        mma_bf16_16816(c[qd], (word << 8) & M2, (word << 10) & M2, (word << 12) & M2,
                       (word << 14) & M2, b[qd].z, b[qd].w);
    }
}

// kModeA: bf16 activations (else int8 from the quantiser).  NT: token
// columns staged (a power of two >= N; columns n >= N repeat token N-1 and
// their results are discarded).
template <bool kModeA, int NT>
__global__ void __launch_bounds__(kThreads, 1)
tl_mma_kernel(const __grid_constant__ GroupArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;                                    // [kWarps][kSlots][2 KB]
    uint4 *xs = reinterpret_cast<uint4 *>(smem + kRingBytes); // staged activations
    __shared__ __align__(8) unsigned long long bars[kWarps][kSlots];
    __shared__ int pend_r[kWarps][kMaxPending];
    __shared__ unsigned long long pend_add[kWarps][kMaxPending];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int v = blockIdx.x * kWarps + warp;
    const int u0 = bnd(a, v), u1 = bnd(a, v + 1);
    const int cu0 = bnd(a, blockIdx.x * kWarps), cu1 = bnd(a, (blockIdx.x + 1) * kWarps);
    const int su = a.R * a.KS;
    const int s_lo = cu0 / su;
    const int n_sl = cu1 > cu0 ? (cu1 - 1) / su - s_lo + 1 : 0;
    const int N = a.N;

    if (threadIdx.x < kWarps * kSlots)
        mbar_init(smem_u32(&bars[0][0]) + 8u * threadIdx.x, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();

    // Weights do not depend on the previous kernel: start the bulk copies
    // before waiting for it.
    const uint32_t ring_w = smem_u32(ring) + warp * (kSlots * kChunkTiles * 512);
    const uint32_t bar_w = smem_u32(&bars[warp][0]);
    Chunk pf;
    pf.seek(a, u0, u1);
    if (lane == 0)
        for (int i = 0; i < kSlots && pf.u < u1; ++i) {
            bulk_load(ring_w + i * (kChunkTiles * 512), pf.src(a), pf.n * 512, bar_w + 8u * i);
            pf.next(a, u1);
        }
    griddep_wait();
    griddep_launch();

    // ---- stage X for this CTA's slices in B-fragment order:
    // word ((((sl*KS + bp)*4 + qd)*NT + n)*4 + t)*4 + w holds x[n'][k], x[n'][k+1],
    // n' = min(n, N-1), k = ((s_lo+sl)*KS + bp)*128 + 16*(2qd + w/2) + 2t + 8*(w%2).
    {
        const int words = n_sl * a.KS * 64 * NT;
        uint32_t *xw = reinterpret_cast<uint32_t *>(xs);
        for (int idx = threadIdx.x; idx < words; idx += kThreads) {
            const int w = idx & 3, tt = (idx >> 2) & 3;
            const int n = min((idx >> 4) % NT, N - 1);
            int rest = (idx >> 4) / NT;
            const int qd = rest & 3;
            rest >>= 2;
            const int bp = rest % a.KS;
            const int sl = rest / a.KS;
            const int k = ((s_lo + sl) * a.KS + bp) * 128 + 16 * (2 * qd + (w >> 1)) + 2 * tt +
                          8 * (w & 1);
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

    // ---- stream the warp's units
    constexpr int XQ = NT * 4;                  // uint4 per 32-column quarter
    constexpr int XB = 4 * XQ;                  // uint4 per 128-column block
    float c[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
    int pend_count = 0;
    int piece_nk = 0;
    Chunk cc;
    cc.seek(a, u0, u1);
    int piece_p = cc.bp == 0 ? 0 : 1;
    int slot = 0;
    uint32_t phases = 0;                        // parity bit per slot
    bool ok = true;

    while (cc.u < u1) {
        const bool got = __all_sync(0xffffffffu, mbar_wait(bar_w + 8u * slot, (phases >> slot) & 1u,
                                                            a.status));
        if (!got) { ok = false; break; }
        phases ^= 1u << slot;
        const uint4 *tiles = reinterpret_cast<const uint4 *>(
            ring + warp * (kSlots * kChunkTiles * 512) + slot * (kChunkTiles * 512)) + lane;
        const uint4 *xb = xs + ((cc.s - s_lo) * a.KS + cc.bp) * XB + (g % NT) * 4 + t;
        if (cc.n == kChunkTiles) {
            // full chunk: load tile i+1 while tile i is multiplied
            uint4 w = tiles[0];
            uint4 b[4];
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) b[qd] = xb[qd * XQ];
#pragma unroll
            for (int i = 0; i < kChunkTiles; ++i) {
                uint4 wn = w, bn[4] = {b[0], b[1], b[2], b[3]};
                if (i + 1 < kChunkTiles) {
                    wn = tiles[(i + 1) * 32];
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd) bn[qd] = xb[(i + 1) * XB + qd * XQ];
                }
                tile_mma(c, w, b);
                w = wn;
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) b[qd] = bn[qd];
            }
        } else {
            for (int i = 0; i < cc.n; ++i) {
                const uint4 w = tiles[i * 32];
                uint4 b[4];
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) b[qd] = xb[i * XB + qd * XQ];
                tile_mma(c, w, b);
            }
        }
        piece_nk += cc.n;
        if (cc.seg_end(a, u1)) {
            // weights decode to +-2: halve (exact)
            pend_count = emit_piece(a, cc.r, cc.s, piece_p, piece_nk, cc.gi, cc.rl, lane,
                                    ((c[0][0] + c[1][0]) + (c[2][0] + c[3][0])) * 0.5f,
                                    ((c[0][1] + c[1][1]) + (c[2][1] + c[3][1])) * 0.5f,
                                    ((c[0][2] + c[1][2]) + (c[2][2] + c[3][2])) * 0.5f,
                                    ((c[0][3] + c[1][3]) + (c[2][3] + c[3][3])) * 0.5f,
                                    pend_r[warp], pend_add[warp], pend_count);
#pragma unroll
            for (int j = 0; j < 4; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
            piece_p = 0;
            piece_nk = 0;
        }
        // refill this slot with the chunk kSlots ahead
        __syncwarp();
        if (lane == 0 && pf.u < u1) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            bulk_load(ring_w + slot * (kChunkTiles * 512), pf.src(a), pf.n * 512, bar_w + 8u * slot);
            pf.next(a, u1);
        }
        cc.next(a, u1);
        slot = slot + 1 == kSlots ? 0 : slot + 1;
    }
    if (!ok) {
        // a copy never landed: drain what is still in flight (bounded), then leave
        for (int i = 0; i < kSlots; ++i) mbar_wait(bar_w + 8u * i, (phases >> i) & 1u, a.status);
        return;
    }
    if (pend_count) commit_pieces(a, pend_r[warp], pend_add[warp], pend_count, lane);
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
                                             (int)(kRingBytes + kSmemLimit)) != cudaSuccess)
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
    int R, KB, KS, S, P;
    long long U, V;
    size_t smem;       // for the given N
    size_t ws_bytes;   // workspace for the given N
};

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// The plan depends on the shapes and the SM count only, never on N, so every
// token is summed in the same order whatever the batch.
void make_plan(const int *Ms, int G, int K, int N, int sms, Plan *p) {
    p->R = 0;
    for (int g = 0; g < G; ++g) p->R += (int)ceil_div(Ms[g], 16);
    p->KB = (int)ceil_div(K, 128);
    p->U = (long long)p->R * p->KB;
    long long ctas = sms;                       // one CTA of kWarps warps per SM
    ctas = std::min<long long>(ctas, ceil_div(p->U, (long long)kWarps * 2));
    if (ctas < 1) ctas = 1;
    p->P = (int)ctas;
    p->V = ctas * kWarps;
    const long long avg = p->U / p->V;
    // Largest slice (in 128-column blocks) that divides KB, keeps every
    // slice segment within two warps (min warp range >= KS - 1) and keeps
    // the staged activations of one CTA within the shared-memory budget at
    // N = 8.  Chosen without looking at N.
    // a CTA covers kWarps consecutive warp ranges of ceil(U/V) units each
    long long cta_units = kWarps * ceil_div(p->U, p->V);
    p->KS = 1;
    for (int d = 1; d <= p->KB && d <= kMaxSlice; ++d) {
        if (p->KB % d != 0 || d > avg + 1) continue;
        const long long su = (long long)p->R * d;
        const long long n_sl = std::min<long long>(p->KB / d, ceil_div(cta_units, su) + 1);
        if ((size_t)n_sl * d * 128 * kNMax * 2 <= kSmemLimit) p->KS = d;
    }
    p->S = p->KB / p->KS;
    if (p->S > kMaxSlices) {                // fewer warps, longer slices
        p->KS = (int)ceil_div(p->KB, kMaxSlices);
        while (p->KB % p->KS) ++p->KS;
        p->S = p->KB / p->KS;
        const long long need_avg = p->KS - 1;       // min warp range >= KS - 1
        long long V = need_avg > 0 ? p->U / need_avg : p->V;
        V = std::max<long long>(kWarps, std::min<long long>(V, p->V)) / kWarps * kWarps;
        p->V = V;
        p->P = (int)(V / kWarps);
    }
    // the per-CTA range may have grown above; size the staging for the final plan
    const long long su = (long long)p->R * p->KS;
    cta_units = kWarps * ceil_div(p->U, p->V);
    const long long n_sl = std::min<long long>(p->S, ceil_div(cta_units, su) + 1);
    const int n = padded_tokens(std::min(std::max(N, 1), kNMax));
    p->smem = (size_t)n_sl * p->KS * 128 * n * 2;
    const size_t cnt_bytes = ((size_t)p->R * 8 + 255) / 256 * 256;
    p->ws_bytes = tl_internal::kStatusBytes + cnt_bytes + (size_t)p->R * p->S * 2 * 16 * n * 4;
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
    make_plan(Ms, G, K, N, sms, &p);
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
    make_plan(Ms, G, K, n, dev.sms, &p);
    if (p.smem > kSmemLimit || p.U >= (1ll << 30)) return TL_ERR_SHAPE;
    if (!ws || ws_bytes < p.ws_bytes) return TL_ERR_WORKSPACE;
    a.R = p.R; a.KB = p.KB; a.KS = p.KS; a.S = p.S; a.K = K; a.U = p.U; a.V = p.V;
    a.L = (int)ceil_div(p.U, p.V);
    const size_t xsz = mode == TL_MODE_BF16 ? 2 : 1;
    a.X = static_cast<const char *>(X) + (size_t)n0 * K * xsz;
    a.s = s ? s + n0 : nullptr;
    a.z = z ? z + n0 : nullptr;
    a.N = n; a.mode = mode; a.out = out;
    const size_t cnt_bytes = ((size_t)p.R * 8 + 255) / 256 * 256;
    char *wsb = static_cast<char *>(ws) + tl_internal::kStatusBytes;
    a.cnt = reinterpret_cast<unsigned long long *>(wsb);
    a.status = static_cast<int *>(ws);
    a.part = reinterpret_cast<float *>(wsb + cnt_bytes);

    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)p.P);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kRingBytes + p.smem;
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
    make_plan(Ms, G, Ws[0].K, kNMax, dev->sms, &p);   // chunks never exceed 8 tokens
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
